"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties one oracle function to an external fact: a published
verification value, a property that characterises linear probing, a library
routine (torch.nn.functional.embedding_bag and its autograd backward,
torch.optim.Adagrad, numpy's float16 cast), a brute-force recomputation, or a
hand-worked example under tests/golden/.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1


# ------------------------------------------------------------------ row-wise Adagrad

def _torch_adagrad(w0, G, acc0, lr, eps):
    p = torch.nn.Parameter(torch.from_numpy(np.asarray(w0, dtype=np.float32).copy()))
    opt = torch.optim.Adagrad([p], lr=lr, eps=eps, initial_accumulator_value=float(acc0))
    p.grad = torch.from_numpy(np.asarray(G, dtype=np.float32))
    opt.step()
    return p.detach().numpy(), opt.state[p]["sum"].numpy()


def test_rowwise_adagrad_one_element_rows_match_torch_adagrad():
    # a row of one element: the row-wise rule is element-wise Adagrad (the library routine)
    rng = np.random.default_rng(31)
    n = 2048
    w0 = rng.uniform(-0.05, 0.05, n).astype(np.float32)
    G = rng.standard_normal(n) * rng.choice([1e-3, 1.0, 30.0], size=n)
    w, acc = oracle.rowwise_adagrad(G, np.arange(n + 1), w0, np.full(n, 0.1, np.float32), 0.01, 1e-8)
    ref_w, ref_acc = _torch_adagrad(w0, G, 0.1, 0.01, 1e-8)
    np.testing.assert_allclose(acc, ref_acc, rtol=2 ** -23, atol=0)
    np.testing.assert_allclose(w, ref_w, rtol=0, atol=2 * np.spacing(np.abs(ref_w)).max())


def test_rowwise_adagrad_equal_gradients_match_elementwise_adagrad():
    # every element of a row with the same gradient g: the row's mean square is g^2, so each
    # element follows torch's element-wise Adagrad from the row's accumulator
    rng = np.random.default_rng(32)
    dims = rng.integers(1, 65, 300)
    goff = np.concatenate([[0], np.cumsum(dims)])
    g_row = rng.standard_normal(dims.size) * 0.5
    G = np.repeat(g_row, dims)
    w0 = rng.uniform(-0.05, 0.05, int(goff[-1])).astype(np.float32)
    w, acc = oracle.rowwise_adagrad(G, goff, w0, np.full(dims.size, 0.1, np.float32), 0.05, 1e-8)
    ref_w, ref_acc = _torch_adagrad(w0, G, 0.1, 0.05, 1e-8)
    # the float32 sum of D equal squares carries up to about D roundings of g^2
    u = 2.0 ** -24
    a_tol = (dims + 2) * u
    np.testing.assert_array_less(np.abs(acc - ref_acc[goff[:-1]]), a_tol * ref_acc[goff[:-1]] + 1e-30)
    step = np.abs(0.05 * G / np.sqrt(np.repeat(ref_acc[goff[:-1]], dims)))
    w_tol = np.repeat(a_tol, dims) * step + 2 * np.spacing(np.abs(ref_w))
    np.testing.assert_array_less(np.abs(w - ref_w), w_tol)


def test_rowwise_adagrad_worked_example_and_order_invariance():
    # hand-worked: g = (1, 7), mean square 25, accumulator 0 -> 25, sqrt 5; lr 5, eps 0:
    # each weight moves by exactly its gradient
    w, acc = oracle.rowwise_adagrad(np.array([1.0, 7.0]), np.array([0, 2]), np.array([10.0, 20.0], np.float32),
                                    np.array([0.0], np.float32), 5.0, 0.0)
    assert np.array_equal(w, np.array([9.0, 13.0], np.float32)) and np.array_equal(acc, np.array([25.0], np.float32))
    # two rows: permuting a row's elements permutes its results (integer gradients: exact sums)
    G = np.array([3.0, -4.0, 12.0, 1.0, 2.0])
    goff = np.array([0, 3, 5])
    w0 = np.array([1.0, 2.0, 3.0, 4.0, 5.0], np.float32)
    a0 = np.array([0.25, 1.5], np.float32)
    w1, a1 = oracle.rowwise_adagrad(G, goff, w0, a0, 0.1, 1e-6)
    perm = np.array([2, 0, 1, 4, 3])
    w2, a2 = oracle.rowwise_adagrad(G[perm], goff, w0[perm], a0, 0.1, 1e-6)
    assert np.array_equal(a1, a2) and np.array_equal(w1[perm], w2)
    assert a1[0] == np.float32(0.25) + np.float32(169.0 / 3) and a1[1] == np.float32(1.5) + np.float32(2.5)
    # half weights: read exactly, rounded to nearest-even like numpy's cast
    wh, _ = oracle.rowwise_adagrad(G, goff, w0.astype(np.float16), a0, 0.1, 1e-6)
    assert np.array_equal(wh, w1.astype(np.float16))


# ------------------------------------------------------------------ fmix64

def _rotl(x, r):
    return ((x << r) | (x >> (64 - r))) & M64


def _murmur3_x64_128(data: bytes, seed: int) -> bytes:
    """MurmurHash3_x64_128 (Appleby), restated from the published algorithm.
    Its finalisation step calls the ORACLE's fmix64, so the verification value
    below pins that function."""
    c1, c2 = 0x87C37B91114253D5, 0x4CF5AD432745937F
    n = len(data)
    h1 = h2 = seed & 0xFFFFFFFF
    nb = n // 16
    for i in range(nb):
        k1 = int.from_bytes(data[16 * i:16 * i + 8], "little")
        k2 = int.from_bytes(data[16 * i + 8:16 * i + 16], "little")
        k1 = (k1 * c1) & M64; k1 = _rotl(k1, 31); k1 = (k1 * c2) & M64; h1 ^= k1
        h1 = _rotl(h1, 27); h1 = (h1 + h2) & M64; h1 = (h1 * 5 + 0x52DCE729) & M64
        k2 = (k2 * c2) & M64; k2 = _rotl(k2, 33); k2 = (k2 * c1) & M64; h2 ^= k2
        h2 = _rotl(h2, 31); h2 = (h2 + h1) & M64; h2 = (h2 * 5 + 0x38495AB5) & M64
    tail = data[16 * nb:]
    k1 = k2 = 0
    for i in range(len(tail) - 1, 7, -1):
        k2 ^= tail[i] << ((i - 8) * 8)
    if len(tail) > 8:
        k2 = (k2 * c2) & M64; k2 = _rotl(k2, 33); k2 = (k2 * c1) & M64; h2 ^= k2
    for i in range(min(len(tail), 8) - 1, -1, -1):
        k1 ^= tail[i] << (i * 8)
    if len(tail) > 0:
        k1 = (k1 * c1) & M64; k1 = _rotl(k1, 31); k1 = (k1 * c2) & M64; h1 ^= k1
    h1 ^= n; h2 ^= n
    h1 = (h1 + h2) & M64; h2 = (h2 + h1) & M64
    h1 = oracle.fmix64(h1); h2 = oracle.fmix64(h2)
    h1 = (h1 + h2) & M64; h2 = (h2 + h1) & M64
    return h1.to_bytes(8, "little") + h2.to_bytes(8, "little")


def test_fmix64_murmur3_verification_value():
    """SMHasher's verification procedure for MurmurHash3_x64_128 yields 0x6384BA69."""
    key = bytes(range(256))
    hashes = b"".join(_murmur3_x64_128(key[:i], 256 - i) for i in range(256))
    final = _murmur3_x64_128(hashes, 0)
    assert int.from_bytes(final[:4], "little") == 0x6384BA69


def test_fmix64_basic_properties():
    assert oracle.fmix64(0) == 0
    rng = np.random.default_rng(1)
    xs = [int(v) for v in rng.integers(0, 2**63, size=2000, dtype=np.int64)]
    assert len({oracle.fmix64(x) for x in xs}) == len(xs)          # injective on a sample
    flips = [bin(oracle.fmix64(x) ^ oracle.fmix64(x ^ 1)).count("1") for x in xs[:500]]
    assert 28 < np.mean(flips) < 36                                  # avalanche


# ------------------------------------------------------------------ table layout

def _tiny_keys(rng, n, n_slots=3):
    raws = rng.choice(1 << 20, size=n, replace=False).astype(np.int64)
    slots = rng.integers(0, n_slots, size=n).astype(np.int64)
    return (slots << 48) | raws


def _home(k, cap):
    return oracle.fmix64(int(k)) & (cap - 1)


@pytest.mark.parametrize("seed,n,cap", [(0, 10, 16), (1, 60, 64), (2, 64, 128), (3, 200, 256), (4, 1, 2)])
def test_layout_characterised_by_linear_probing(seed, n, cap):
    """Every key sits at the first slot of its cyclic probe path that no EARLIER
    key took: all slots between its home and its slot hold earlier keys."""
    rng = np.random.default_rng(seed)
    keys = _tiny_keys(rng, n)
    T = oracle.Table(keys, cap, [4, 4, 4])
    sk, sr = T.layout()
    pos = {int(k): i for i, k in enumerate(keys)}
    occupied = np.nonzero(sk != -1)[0]
    assert len(occupied) == n and sorted(sk[occupied].tolist()) == sorted(keys.tolist())
    max_probe = 0
    for p in occupied:
        k = int(sk[p])
        assert sr[p] == pos[k]
        h = _home(k, cap)
        d = (p - h) % cap
        for j in range(d):
            q = (h + j) % cap
            assert sk[q] != -1 and pos[int(sk[q])] < pos[k]
        max_probe = max(max_probe, d + 1)
    assert T.max_probe == max_probe
    # longest cyclic run of occupied slots, counted directly
    occ = np.concatenate([sk != -1, sk != -1])
    best = run = 0
    for o in occ:
        run = run + 1 if o else 0
        best = max(best, run)
    assert T.max_cluster == min(best, cap)


def test_layout_occupied_set_independent_of_insert_order():
    rng = np.random.default_rng(7)
    keys = _tiny_keys(rng, 500)
    a, _ = oracle.Table(keys, 1024, [4, 4, 4]).layout()
    b, _ = oracle.Table(keys[rng.permutation(500)], 1024, [4, 4, 4]).layout()
    assert np.array_equal(a != -1, b != -1)
    assert not np.array_equal(a, b)    # assignment does depend on the order


def test_resolve_brute_force():
    rng = np.random.default_rng(3)
    keys = _tiny_keys(rng, 100)
    T = oracle.Table(keys, 256, [4, 4, 4])
    sk, _ = T.layout()
    absent = _tiny_keys(np.random.default_rng(99), 200)
    absent = absent[~np.isin(absent, keys)]
    q = np.concatenate([keys, absent, [-1]])
    slot, row = T.resolve(q)
    for i, k in enumerate(q):
        where = np.nonzero(sk == k)[0] if k != -1 else []
        if len(where):
            assert slot[i] == where[0] and keys[row[i]] == k
        else:
            assert slot[i] == -1 and row[i] == -1


def test_build_rejects_bad_tables():
    with pytest.raises(oracle.OracleError, match="duplicate"):
        oracle.Table(np.array([1, 2, 1]), 8, [4])
    with pytest.raises(oracle.OracleError, match="reserved"):
        oracle.Table(np.array([1, -1]), 8, [4])
    with pytest.raises(oracle.OracleError, match="bad slot"):
        oracle.Table(np.array([(3 << 48) | 1]), 8, [4, 4])
    with pytest.raises(oracle.OracleError, match="invalid"):
        oracle.Table(np.array([1, 2]), 6, [4])


# ------------------------------------------------------------------ golden fixtures

def test_golden_key_layout():
    g = json.load(open(os.path.join(GOLDEN, "unified_key_layout.json")))
    for c in g["cases"]:
        k = c["key"]
        assert (c["slot"] << 48) | c["raw"] == k
        # the oracle reads the slot field from the high 16 bits: a table whose
        # slots have distinct dims places the row accordingly
        dims = [1] * 32768
        dims[c["slot"]] = 3
        T = oracle.Table(np.array([k], dtype=np.int64), 2, dims)
        assert T.elem_offsets().tolist() == [0, 3]


def test_golden_csr_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "csr_worked_example.json")))
    T = oracle.Table(np.array(g["table_keys"], dtype=np.int64), g["capacity"], g["dims"])
    values = np.array(g["values"], dtype=np.float32).reshape(-1)
    off = np.array(g["offsets"]); keys = np.array(g["keys"], dtype=np.int64)
    grad = np.array(g["grad_out"], dtype=np.float32)
    for pool in ("sum", "mean"):
        out, _ = T.forward(off, keys, pool, "f32", values)
        np.testing.assert_allclose(out, np.array(g[pool]), rtol=1e-15, atol=0)
        uk, _, goff, G, _ = T.backward(off, keys, pool, grad)
        assert uk.tolist() == g["unique_keys"]
        for i, k in enumerate(uk):
            np.testing.assert_allclose(G[goff[i]:goff[i + 1]], g["G_" + pool][str(int(k))], rtol=1e-15)


# ------------------------------------------------------------------ pooling vs torch EmbeddingBag

def _random_case(seed, n_keys=300, n_slots=3, D=8, B=40, max_len=12, absent_p=0.2, wd=np.float32):
    rng = np.random.default_rng(seed)
    keys = np.empty(0, dtype=np.int64)
    per = n_keys // n_slots
    for s in range(n_slots):
        keys = np.concatenate([keys, (np.int64(s) << 48) | rng.choice(1 << 30, size=per, replace=False)])
    keys = keys[rng.permutation(keys.size)]
    values = rng.standard_normal((keys.size, D)).astype(wd)
    L = rng.integers(0, max_len + 1, size=B * n_slots)
    off = np.concatenate([[0], np.cumsum(L)])
    q = np.empty(off[-1], dtype=np.int64)
    for bag in range(B * n_slots):
        s = bag % n_slots
        mine = keys[(keys >> 48) == s]
        pick = mine[rng.integers(0, mine.size, size=L[bag])]
        miss = rng.random(L[bag]) < absent_p
        pick[miss] = (np.int64(s) << 48) | ((1 << 31) + rng.integers(0, 1000, size=miss.sum()))
        q[off[bag]:off[bag + 1]] = pick
    grad = rng.standard_normal((B, n_slots * D)).astype(np.float32)
    return keys, values, off, q, grad


@pytest.mark.parametrize("wd", [np.float32, np.float16], ids=["f32", "f16"])
@pytest.mark.parametrize("pool", ["sum", "mean"])
def test_forward_matches_torch_embedding_bag(pool, wd):
    """Float32 and float16 rows: the half rows are read by the oracle's own
    half loader and by numpy's exact half -> double conversion here, so a
    wrong element width, offset or conversion in the former fails."""
    keys, values, off, q, _ = _random_case(11, absent_p=0.0, wd=wd)
    n_slots, D = 3, 8
    T = oracle.Table(keys, 1024, [D] * n_slots)
    out, A = T.forward(off, q, pool, "f16" if wd == np.float16 else "f32", values.reshape(-1))
    # library routine: EmbeddingBag over dense row indices (independent dict lookup)
    idx = {int(k): i for i, k in enumerate(keys)}
    flat = torch.tensor([idx[int(k)] for k in q], dtype=torch.int64)
    ref = torch.nn.functional.embedding_bag(flat, torch.from_numpy(values.astype(np.float64)),
                                            torch.from_numpy(off[:-1]), mode=pool)
    np.testing.assert_allclose(out.reshape(-1, D), ref.numpy(), rtol=1e-13, atol=1e-13)
    assert np.all(A.reshape(-1, D) >= np.abs(out.reshape(-1, D)) - 1e-12)


@pytest.mark.parametrize("pool", ["sum", "mean"])
def test_backward_matches_torch_autograd(pool):
    keys, values, off, q, grad = _random_case(12, absent_p=0.0)
    n_slots, D = 3, 8
    T = oracle.Table(keys, 1024, [D] * n_slots)
    uk, rows, goff, G, _ = T.backward(off, q, pool, grad)
    idx = {int(k): i for i, k in enumerate(keys)}
    flat = torch.tensor([idx[int(k)] for k in q], dtype=torch.int64)
    W = torch.from_numpy(values).double().requires_grad_(True)
    y = torch.nn.functional.embedding_bag(flat, W, torch.from_numpy(off[:-1]), mode=pool)
    # pooled rows are bags in sample-major order: bag b*S+s <- grad_out[b, s*D:(s+1)*D]
    y.backward(torch.from_numpy(grad).double().reshape(-1, D))
    ref = W.grad.numpy()
    assert set(uk.tolist()) == set(q.tolist())
    assert sorted(rows.tolist()) == sorted(np.nonzero(np.abs(ref).sum(1) > 0)[0].tolist())
    for i, r in enumerate(rows):
        np.testing.assert_allclose(G[goff[i]:goff[i + 1]], ref[r], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("wd", [np.float32, np.float16], ids=["f32", "f16"])
def test_pooling_brute_force_with_misses_and_special_cases(wd):
    keys, values, off, q, grad = _random_case(13, absent_p=0.3, max_len=6, wd=wd)
    n_slots, D = 3, 8
    T = oracle.Table(keys, 1024, [D] * n_slots)
    table = {int(k): values[i].astype(np.float64) for i, k in enumerate(keys)}
    wname = "f16" if wd == np.float16 else "f32"
    s_out, _ = T.forward(off, q, "sum", wname, values.reshape(-1))
    m_out, _ = T.forward(off, q, "mean", wname, values.reshape(-1))
    s_out = s_out.reshape(-1, D); m_out = m_out.reshape(-1, D)
    for bag in range(off.size - 1):
        ks = q[off[bag]:off[bag + 1]]
        hits = [table[int(k)] for k in ks if int(k) in table]
        exp = np.array([math.fsum(h[j] for h in hits) for j in range(D)]) if hits else np.zeros(D)
        np.testing.assert_allclose(s_out[bag], exp, rtol=1e-13, atol=1e-13)
        L = ks.size
        if L == 0 or not hits:
            assert np.all(s_out[bag] == 0) and np.all(m_out[bag] == 0)      # all-miss / empty bag -> 0
        else:
            np.testing.assert_array_equal(m_out[bag], s_out[bag] / L)        # mean == sum / L
        if L == 1 and hits:
            np.testing.assert_array_equal(s_out[bag], hits[0])               # L=1 sum is the row


def test_backward_brute_force_and_single_hit():
    keys, values, off, q, grad = _random_case(14, absent_p=0.25)
    n_slots, D = 3, 8
    T = oracle.Table(keys, 1024, [D] * n_slots)
    present = set(int(k) for k in keys)
    for pool in ("sum", "mean"):
        uk, rows, goff, G, A = T.backward(off, q, pool, grad)
        contrib = {}
        for bag in range(off.size - 1):
            L = off[bag + 1] - off[bag]
            for k in q[off[bag]:off[bag + 1]]:
                if int(k) in present:
                    b, s = divmod(bag, n_slots)
                    contrib.setdefault(int(k), []).append(
                        grad[b, s * D:(s + 1) * D].astype(np.float64) * (1.0 / L if pool == "mean" else 1.0))
        assert uk.tolist() == sorted(contrib)
        for i, k in enumerate(uk):
            terms = contrib[int(k)]
            exp = [math.fsum(t[j] for t in terms) for j in range(D)]
            np.testing.assert_allclose(G[goff[i]:goff[i + 1]], exp, rtol=1e-13, atol=1e-13)
            if len(terms) == 1:
                np.testing.assert_array_equal(G[goff[i]:goff[i + 1]], terms[0])
            np.testing.assert_allclose(A[goff[i]:goff[i + 1]],
                                       [math.fsum(abs(t[j]) for t in terms) for j in range(D)], rtol=1e-13)


def test_ragged_dims_offsets_and_pooling():
    rng = np.random.default_rng(5)
    dims = [8, 16, 4]
    keys = np.concatenate([(np.int64(s) << 48) | rng.choice(1 << 20, size=20, replace=False) for s in range(3)])
    keys = keys[rng.permutation(keys.size)]
    T = oracle.Table(keys, 128, dims)
    off_e = T.elem_offsets()
    d = np.array([dims[k >> 48] for k in keys])
    assert off_e.tolist() == [0] + np.cumsum(d).tolist()
    values = rng.standard_normal(off_e[-1]).astype(np.float32)
    # one sample, one bag per slot, each bag pooling every key of its slot
    bags = [keys[(keys >> 48) == s] for s in range(3)]
    off = np.array([0] + np.cumsum([b.size for b in bags]).tolist())
    out, _ = T.forward(off, np.concatenate(bags), "sum", "f32", values)
    pos = {int(k): i for i, k in enumerate(keys)}
    exp = np.concatenate([
        np.sum([values[off_e[pos[int(k)]]:off_e[pos[int(k)] + 1]].astype(np.float64) for k in bags[s]], axis=0)
        for s in range(3)])
    np.testing.assert_allclose(out.reshape(-1), exp, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ Adagrad

@pytest.mark.parametrize("wd", [np.float32, np.float16])
def test_adagrad_matches_torch_optim_adagrad(wd):
    rng = np.random.default_rng(21)
    n = 4096
    w0 = (rng.uniform(-0.05, 0.05, n)).astype(wd)
    acc0 = np.full(n, 0.1, dtype=np.float32)
    G = rng.standard_normal(n) * rng.choice([1e-3, 1.0, 30.0], size=n)
    G[:64] = 0.0
    lr, eps = 0.01, 1e-8
    w, acc = oracle.adagrad(G, w0, acc0, lr, eps)
    # library routine: torch.optim.Adagrad, float32, initial accumulator 0.1
    p = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float32)))
    opt = torch.optim.Adagrad([p], lr=lr, eps=eps, initial_accumulator_value=0.1)
    p.grad = torch.from_numpy(G.astype(np.float32))
    opt.step()
    ref_w = p.detach().numpy().astype(wd)
    ref_acc = opt.state[p]["sum"].numpy()
    np.testing.assert_allclose(acc, ref_acc, rtol=2 ** -23, atol=0)
    if wd == np.float32:
        np.testing.assert_allclose(w, ref_w, rtol=0, atol=2 * np.spacing(np.abs(ref_w)).max())
    else:
        # half results may differ only where float32 noise straddles a rounding boundary
        assert np.mean(w == ref_w) > 0.999
        np.testing.assert_allclose(w.astype(np.float32), ref_w.astype(np.float32), rtol=0,
                                   atol=float(np.spacing(np.float16(0.06))))
    # g = 0 leaves the row bit-identical (features absent from a batch are untouched)
    assert np.array_equal(w[:64], w0[:64]) and np.array_equal(acc[:64], acc0[:64])


def test_adagrad_single_hit_closed_form():
    rng = np.random.default_rng(22)
    n = 2000
    w0 = rng.uniform(-0.05, 0.05, n).astype(np.float32)
    acc0 = rng.uniform(0.01, 2.0, n).astype(np.float32)
    g = rng.standard_normal(n).astype(np.float32).astype(np.float64)
    lr, eps = 0.01, 1e-8
    w, acc = oracle.adagrad(g, w0, acc0, lr, eps)
    acc_cf = acc0.astype(np.float64) + g * g
    w_cf = w0.astype(np.float64) - lr * g / (np.sqrt(acc_cf) + eps)
    np.testing.assert_allclose(acc, acc_cf, rtol=3e-7)
    np.testing.assert_allclose(w, w_cf, rtol=0, atol=4 * np.spacing(np.float32(0.06)))


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(23)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 0.05,
        rng.standard_normal(2000).astype(np.float32) * 1e-6,          # subnormal halves
        np.float32([65504, 65520, 65519.99, 1e9, -1e9, 0.0, -0.0, 6e-8, 3e-8, np.inf, -np.inf]),
    ])
    # exact halfway cases between adjacent halves
    h = rng.integers(0, 0x7BFF, size=2000, dtype=np.uint16).view(np.float16)
    mid = ((h.astype(np.float64) + np.nextafter(h, np.float16(np.inf)).astype(np.float64)) / 2).astype(np.float32)
    x = np.concatenate([x, mid])
    assert np.array_equal(oracle.f32_to_f16_bits(x), x.astype(np.float16).view(np.uint16))


def test_master_copy_rows_are_the_masters_rounded_to_nearest_even():
    rng = np.random.default_rng(7)
    m = np.concatenate([rng.uniform(-0.05, 0.05, 4096).astype(np.float32),
                        # exact ties between neighbouring halves go to the even one
                        np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, -(1 + 2.0 ** -11), 65504.0, 1e-8],
                                 dtype=np.float32)])
    c = oracle.f16_copy(m)
    assert c.dtype == np.float16
    assert np.array_equal(c.view(np.uint16), m.astype(np.float16).view(np.uint16))
    assert c[-5] == np.float16(1.0) and c[-4] == np.float16(1 + 2.0 ** -9) and c[-3] == np.float16(-1.0)



# ------------------------------------------------------------------ FTRL-Proximal

def test_ftrl_without_regularisation_is_adagrad():
    """With lambda1 = lambda2 = 0, FTRL-Proximal with per-coordinate rates
    eta_t = alpha / (beta + sqrt(n_t)) is online gradient descent with those
    rates (McMahan et al., KDD 2013, section 3.1: the FTRL-Proximal and OGD
    updates coincide), i.e. Adagrad with lr = alpha and eps = beta, provided
    the starting weight is the one z encodes, w_0 = -eta_0 z_0.  So several
    oracle FTRL steps must follow torch.optim.Adagrad (float64) from that start.
    A wrong sign, a dropped sigma * w term, or sqrt(n) taken before instead of
    after the update breaks the agreement."""
    rng = np.random.default_rng(21)
    m, alpha, beta, n0 = 4000, 0.05, 0.7, 0.1
    w0 = rng.uniform(-0.05, 0.05, m).astype(np.float32)
    z = (-w0.astype(np.float64) * (beta + math.sqrt(n0)) / alpha).astype(np.float32)
    n = np.full(m, n0, np.float32)
    w = w0.copy()
    p = torch.from_numpy(w0.astype(np.float64)).requires_grad_(True)
    opt = torch.optim.Adagrad([p], lr=alpha, eps=beta, initial_accumulator_value=n0)
    for step in range(6):
        g = rng.standard_normal(m) * (0.3 if step % 2 else 2.0)
        w, n, z = oracle.ftrl(g, w, n, z, alpha, beta, 0.0, 0.0)
        p.grad = torch.from_numpy(g.astype(np.float32).astype(np.float64))
        opt.step()
        ref = p.detach().numpy()
        np.testing.assert_allclose(w, ref, rtol=2e-5, atol=2e-5 * np.abs(ref).max())


def test_ftrl_weight_is_the_proximal_minimiser():
    """The closed-form weight is the minimiser of the per-coordinate objective
    z w + lambda1 |w| + (1/2) ((beta + sqrt(n)) / alpha + lambda2) w^2
    (McMahan et al. 2013, Algorithm 1 and its derivation); checked against a
    numerical minimisation, which pins the signs and where lambda1 and
    lambda2 enter.  One step from w = 0 (so z' = z + g exactly)."""
    from scipy.optimize import minimize_scalar
    rng = np.random.default_rng(22)
    alpha, beta, l1, l2 = 0.1, 1.0, 0.4, 0.3
    m = 300
    g = rng.standard_normal(m) * 1.5
    w, n, z = oracle.ftrl(g, np.zeros(m, np.float32), np.full(m, 0.25, np.float32),
                          rng.standard_normal(m).astype(np.float32), alpha, beta, l1, l2)
    zeros = 0
    for i in range(m):
        q = (beta + math.sqrt(float(n[i]))) / alpha + l2
        f = lambda x: float(z[i]) * x + l1 * abs(x) + 0.5 * q * x * x
        r = minimize_scalar(f, bounds=(-50.0, 50.0), method="bounded", options={"xatol": 1e-12})
        assert abs(float(w[i]) - r.x) <= 1e-6 * max(1.0, abs(r.x)), (i, w[i], r.x)
        zeros += w[i] == 0
    assert 0 < zeros < m                         # both branches exercised


def test_ftrl_state_invariants():
    """n accumulates g^2 exactly as the Adagrad accumulator does (same float32
    operations); with w = 0 the z update is z + g; lambda1 above every |z|
    makes every weight exactly 0 (the sparsity FTRL-Proximal is used for)."""
    rng = np.random.default_rng(23)
    m = 1000
    G = rng.standard_normal(m)
    w0 = rng.uniform(-0.05, 0.05, m).astype(np.float32)
    n0 = np.full(m, 0.1, np.float32)
    z0 = rng.standard_normal(m).astype(np.float32)
    _, n1, _ = oracle.ftrl(G, w0, n0, z0, 0.05, 1.0, 0.0, 0.0)
    _, acc1 = oracle.adagrad(G, w0, n0, 0.05, 1e-8)
    assert np.array_equal(n1.view(np.uint32), acc1.view(np.uint32))
    _, _, z1 = oracle.ftrl(G, np.zeros(m, np.float32), n0, z0, 0.05, 1.0, 0.0, 0.0)
    assert np.array_equal(z1, (z0 + G.astype(np.float32)).astype(np.float32))
    wbig, _, _ = oracle.ftrl(G, w0, n0, z0, 0.05, 1.0, 1e6, 0.0)
    assert np.all(wbig == 0)
    wh, _, _ = oracle.ftrl(G, w0.astype(np.float16), n0, z0, 0.05, 1.0, 0.1, 0.2)
    wf, _, _ = oracle.ftrl(G, w0.astype(np.float16).astype(np.float32), n0, z0, 0.05, 1.0, 0.1, 0.2)
    assert wh.dtype == np.float16 and np.array_equal(wh, wf.astype(np.float16))   # half: read exactly, RNE out
