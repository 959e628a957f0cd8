"""Seeded synthetic inputs for the unified-hash-table embedding step.

Input generation only: this module builds keys, CSR batches, initial weights,
initial accumulators and upstream gradients.  It holds none of the step's own
arithmetic (no hashing of keys into the table, no probing, no pooling, no
gradient reduction, no optimizer); both the CUDA path and the oracle consume
the arrays it returns.

Every random number is a pure function of (seed, stream, counter): a
splitmix64-style mixer (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014, the SplitMix64 output function) applied to a
64-bit counter.  It is written with wrapping int64 torch ops, so the same call
gives the same integers on the CPU and on a CUDA device.  Draws that go through
transcendental functions (the Box-Muller normals for ``grad_out``) may differ
in the last bit between devices; parity always feeds ONE generated array to
both sides, so that never matters.

Workload recipe (the five configurations of the embedding-step benchmark):

* keys: ``key = (slot << 48) | raw`` (unified hash table key layout: low 48
  bits raw feature id, high 16 bits table id; Tencent PCG DataFun talk,
  "计算优化" paragraph on the Unified Hash Table).  Per slot ``s`` the table
  holds ranks ``0..V_s-1``; ``raw = (a_s * rank + c_s) mod 2^48`` with an odd
  seeded ``a_s`` (a bijection, so raws never collide).
* keys-array order (the order handed to table creation) is a seeded
  pseudo-random permutation of all (slot, rank) pairs, so hot rows carry no
  artificial locality.
* bags: ``B * S`` bags in sample-major order (bag = b * S + s).  Lengths from
  the configuration's distribution; ids Zipf(s) over ranks of the bag's slot
  (weight ``(rank + 1) ** -s``), drawn by inverse CDF on a float64 table.
* absent keys: with probability ``absent`` an occurrence takes rank
  ``V_s + rank`` instead, which is never in the table (same Zipf popularity).
* initial weights ``U(-0.05, 0.05)`` per element (float32, then float16 for
  half tables); initial accumulators the constant ``acc0``; ``grad_out``
  ``N(0, grad_std^2)`` per element, float32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

__all__ = [
    "Config", "CONFIGS", "config", "scaled",
    "mix64", "uniform01",
    "table_keys", "batch", "w0_values", "w0_rows", "grad_out", "elem_offsets",
    "Workload", "make",
]

_M64 = (1 << 64) - 1


def _s64(c: int) -> int:
    """An unsigned 64-bit constant as the signed int64 torch stores."""
    c &= _M64
    return c - (1 << 64) if c >= (1 << 63) else c


_GOLDEN = _s64(0x9E3779B97F4A7C15)
_MUL1 = _s64(0xBF58476D1CE4E5B9)
_MUL2 = _s64(0x94D049BB133111EB)
_SEEDMUL = _s64(0xD1B54A32D192ED03)
_STREAMMUL = _s64(0xAEF17502108EF2D9)

# purpose streams: one independent sub-stream per kind of draw
STREAM = {
    "vocab": 1, "affine": 2, "order": 3, "len": 4, "id": 5, "absent": 6,
    "w0": 7, "g1": 8, "g2": 9,
}


def _lsr(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def mix64(seed: int, stream: int, counter: torch.Tensor) -> torch.Tensor:
    """SplitMix64 output function of ``seed*A + stream*B + counter`` (wrapping)."""
    x = counter.to(torch.int64) + _s64(seed * _SEEDMUL + stream * _STREAMMUL + _GOLDEN)
    x = (x ^ _lsr(x, 30)) * _MUL1
    x = (x ^ _lsr(x, 27)) * _MUL2
    return x ^ _lsr(x, 31)


def uniform01(seed: int, stream: int, counter: torch.Tensor) -> torch.Tensor:
    """float64 in [0, 1): the top 53 bits of the mixed counter."""
    return _lsr(mix64(seed, stream, counter), 11).to(torch.float64) * (2.0 ** -53)


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    n_slots: int
    vocab: Tuple[int, ...]          # keys per slot, V_s
    dims: Tuple[int, ...]           # embedding dim per slot
    wdtype: str                     # "f32" | "f16" | "f16m" (f32 master + f16 copy; accumulator always f32)
    batch: int                      # samples B; bags = B * n_slots
    bag_len: Tuple                  # ("uniform", lo, hi) | ("geometric", p, cap) | ("zipf", s, lo, hi)
    zipf_s: float
    absent: float
    pool: str                       # "sum" | "mean"
    lr: float
    eps: float
    acc0: float
    grad_std: float
    seed: int = 0

    @property
    def n_keys(self) -> int:
        return int(sum(self.vocab))

    @property
    def n_bags(self) -> int:
        return self.batch * self.n_slots

    @property
    def sum_dims(self) -> int:
        return int(sum(self.dims))

    @property
    def capacity(self) -> int:
        """Smallest power of two holding the keys at load factor <= 0.5."""
        c = 1
        while c < 2 * self.n_keys:
            c <<= 1
        return c

    @property
    def uniform_dim(self) -> bool:
        return len(set(self.dims)) == 1


def _log_uniform_vocab(seed: int, n_slots: int, lo: float, hi: float, total: int) -> Tuple[int, ...]:
    u = uniform01(seed, STREAM["vocab"], torch.arange(n_slots)).numpy()
    v = np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    v = np.rint(v * (total / v.sum())).astype(np.int64)
    v[-1] += total - int(v.sum())
    return tuple(int(x) for x in v)


def _make_configs() -> Dict[int, Config]:
    c = {}
    c[1] = Config("tiny-4slot-16d-f32", 4, (16384,) * 4, (16,) * 4, "f32", 256,
                  ("uniform", 1, 8), 1.05, 0.0, "sum", 0.01, 1e-8, 0.1, 1.0)
    c[2] = Config("26slot-10M-64d-f32-mean", 26, _log_uniform_vocab(0, 26, 1e3, 2e6, 10_000_000),
                  (64,) * 26, "f32", 16384, ("uniform", 1, 20), 1.1, 0.02, "mean", 0.05, 1e-8, 0.1, 1.0)
    c[3] = Config("100slot-50M-32d-f16", 100, (500_000,) * 100, (32,) * 100, "f16", 65536,
                  ("uniform", 1, 10), 1.2, 0.0, "sum", 0.01, 1e-6, 0.1, 1.0)
    c[4] = Config("40slot-20M-ragged-f32", 40, (500_000,) * 40,
                  tuple((8, 16, 32, 64, 128)[s % 5] for s in range(40)), "f32", 32768,
                  ("geometric", 0.2, 64), 1.05, 0.0, "sum", 0.02, 1e-8, 0.1, 1.0)
    c[5] = Config("large-64slot-100M-128d-f16-mean", 64, (1_562_500,) * 64, (128,) * 64, "f16", 131072,
                  ("zipf", 1.1, 1, 256), 1.1, 0.05, "mean", 0.01, 1e-8, 0.1, 0.1)
    return c


CONFIGS: Dict[int, Config] = _make_configs()


def config(i: int) -> Config:
    return CONFIGS[i]


def scaled(cfg: Config, vocab_div: int = 1, batch_div: int = 1, name: Optional[str] = None,
           **override) -> Config:
    """A smaller copy of a configuration with the same structure."""
    vocab = tuple(max(8, v // vocab_div) for v in cfg.vocab)
    fields = dict(vocab=vocab, batch=max(1, cfg.batch // batch_div),
                  name=name or f"{cfg.name}/v{vocab_div}b{batch_div}")
    fields.update(override)
    return dataclasses.replace(cfg, **fields)


# ---------------------------------------------------------------- keys

def _slot_affine(cfg: Config, dev) -> Tuple[torch.Tensor, torch.Tensor]:
    s = torch.arange(cfg.n_slots, device=dev)
    a = (_lsr(mix64(cfg.seed, STREAM["affine"], 2 * s), 16)) | 1          # odd, < 2^48
    c = _lsr(mix64(cfg.seed, STREAM["affine"], 2 * s + 1), 16)             # < 2^48
    return a, c


def _raw(a: torch.Tensor, c: torch.Tensor, rank: torch.Tensor) -> torch.Tensor:
    return (a * rank + c) & ((1 << 48) - 1)


def table_keys(cfg: Config, device="cpu") -> torch.Tensor:
    """int64[N] keys in keys-array order (the order given to table creation)."""
    dev = torch.device(device)
    V = torch.tensor(cfg.vocab, dtype=torch.int64, device=dev)
    base = torch.cumsum(V, 0) - V
    n = cfg.n_keys
    gid = torch.arange(n, dtype=torch.int64, device=dev)
    slot = torch.repeat_interleave(torch.arange(cfg.n_slots, device=dev), V)
    rank = gid - base[slot]
    a, c = _slot_affine(cfg, dev)
    keys = (slot << 48) | _raw(a[slot], c[slot], rank)
    del rank, gid
    # seeded permutation: sort by a bijective hash of the global index (no ties)
    order = torch.argsort(mix64(cfg.seed, STREAM["order"], torch.arange(n, device=dev)))
    return keys[order].contiguous()


# ---------------------------------------------------------------- batches

def _len_cdf(cfg: Config) -> Tuple[np.ndarray, int]:
    kind = cfg.bag_len[0]
    if kind == "geometric":
        p, cap = cfg.bag_len[1], cfg.bag_len[2]
        k = np.arange(1, cap + 1, dtype=np.float64)
        pmf = (1.0 - p) ** (k - 1) * p
        cdf = np.cumsum(pmf)
        cdf[-1] = np.inf  # the cap absorbs the tail
        return cdf, 1
    if kind == "zipf":
        s, lo, hi = cfg.bag_len[1], cfg.bag_len[2], cfg.bag_len[3]
        k = np.arange(lo, hi + 1, dtype=np.float64)
        w = k ** -s
        cdf = np.cumsum(w) / w.sum()
        cdf[-1] = np.inf
        return cdf, lo
    raise ValueError(kind)


def _zipf_cdf(V: int, s: float) -> np.ndarray:
    w = np.arange(1, V + 1, dtype=np.float64) ** -s
    cdf = np.cumsum(w) / w.sum()
    cdf[-1] = np.inf
    return cdf


def bag_lengths(cfg: Config, device="cpu") -> torch.Tensor:
    dev = torch.device(device)
    q = torch.arange(cfg.n_bags, dtype=torch.int64, device=dev)
    u = uniform01(cfg.seed, STREAM["len"], q)
    if cfg.bag_len[0] == "uniform":
        lo, hi = cfg.bag_len[1], cfg.bag_len[2]
        return lo + torch.floor(u * (hi - lo + 1)).to(torch.int64)
    cdf, lo = _len_cdf(cfg)
    return lo + torch.searchsorted(torch.from_numpy(cdf).to(dev), u, right=True)


def batch(cfg: Config, device="cpu") -> Tuple[torch.Tensor, torch.Tensor]:
    """(offsets int64[B*S+1], keys int64[nnz]) in CSR, bag = b * S + s."""
    dev = torch.device(device)
    L = bag_lengths(cfg, dev)
    offsets = torch.zeros(cfg.n_bags + 1, dtype=torch.int64, device=dev)
    torch.cumsum(L, 0, out=offsets[1:])
    nnz = int(offsets[-1])
    slot = torch.repeat_interleave(torch.arange(cfg.n_bags, device=dev) % cfg.n_slots, L)
    del L
    occ = torch.arange(nnz, dtype=torch.int64, device=dev)
    u = uniform01(cfg.seed, STREAM["id"], occ)
    rank = torch.empty(nnz, dtype=torch.int64, device=dev)
    by_v: Dict[int, List[int]] = {}
    for s, v in enumerate(cfg.vocab):
        by_v.setdefault(v, []).append(s)
    for v, slots in by_v.items():
        cdf = torch.from_numpy(_zipf_cdf(v, cfg.zipf_s)).to(dev)
        if len(by_v) == 1:
            rank = torch.searchsorted(cdf, u, right=True)
        else:
            m = torch.isin(slot, torch.tensor(slots, device=dev))
            rank[m] = torch.searchsorted(cdf, u[m], right=True)
    del u
    if cfg.absent > 0:
        ua = uniform01(cfg.seed, STREAM["absent"], occ)
        V = torch.tensor(cfg.vocab, dtype=torch.int64, device=dev)
        rank = torch.where(ua < cfg.absent, rank + V[slot], rank)
        del ua
    a, c = _slot_affine(cfg, dev)
    keys = (slot << 48) | _raw(a[slot], c[slot], rank)
    return offsets, keys.contiguous()


# ---------------------------------------------------------------- values

def elem_offsets(cfg: Config, keys: torch.Tensor) -> torch.Tensor:
    """int64[N+1] element offset of each keys-array row in the ragged values array."""
    dims = torch.tensor(cfg.dims, dtype=torch.int64, device=keys.device)
    d = dims[keys >> 48]
    off = torch.zeros(keys.numel() + 1, dtype=torch.int64, device=keys.device)
    torch.cumsum(d, 0, out=off[1:])
    return off


def _w0_from_elem(cfg: Config, e: torch.Tensor) -> torch.Tensor:
    w = (-0.05 + 0.1 * uniform01(cfg.seed, STREAM["w0"], e)).to(torch.float32)
    return w.to(torch.float16) if cfg.wdtype == "f16" else w


def w0_values(cfg: Config, n_elems: int, device="cpu", chunk: int = 1 << 28,
              out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Initial weights for the whole ragged values array (keys-array row order)."""
    dev = torch.device(device)
    dt = torch.float16 if cfg.wdtype == "f16" else torch.float32
    if out is None:
        out = torch.empty(n_elems, dtype=dt, device=dev)
    for s in range(0, n_elems, chunk):
        e = torch.arange(s, min(n_elems, s + chunk), dtype=torch.int64, device=dev)
        out[s:s + e.numel()] = _w0_from_elem(cfg, e)
    return out


def w0_rows(cfg: Config, elem_off: torch.Tensor, rows: torch.Tensor, dims_of_rows: torch.Tensor):
    """Initial weights of selected keys-array rows, concatenated (ragged)."""
    if rows.numel() == 0:
        return _w0_from_elem(cfg, torch.zeros(0, dtype=torch.int64))
    start = elem_off[rows]
    rep = torch.repeat_interleave(start, dims_of_rows)
    within = torch.arange(int(dims_of_rows.sum()), dtype=torch.int64) - \
        torch.repeat_interleave(torch.cumsum(dims_of_rows, 0) - dims_of_rows, dims_of_rows)
    return _w0_from_elem(cfg, rep + within)


def grad_out(cfg: Config, device="cpu", chunk: int = 1 << 27) -> torch.Tensor:
    """float32[B, sum(dims)] upstream gradient of the pooled output."""
    dev = torch.device(device)
    n = cfg.batch * cfg.sum_dims
    out = torch.empty(n, dtype=torch.float32, device=dev)
    for s in range(0, n, chunk):
        e = torch.arange(s, min(n, s + chunk), dtype=torch.int64, device=dev)
        u1 = uniform01(cfg.seed, STREAM["g1"], e)
        u2 = uniform01(cfg.seed, STREAM["g2"], e)
        z = torch.sqrt(-2.0 * torch.log1p(-u1)) * torch.cos((2.0 * math.pi) * u2)
        out[s:s + e.numel()] = (cfg.grad_std * z).to(torch.float32)
    return out.view(cfg.batch, cfg.sum_dims)


@dataclasses.dataclass
class Workload:
    cfg: Config
    keys: torch.Tensor          # table keys, keys-array order
    offsets: torch.Tensor       # CSR offsets over bags
    qkeys: torch.Tensor         # CSR keys (occurrences)
    values: Optional[torch.Tensor]
    grad: torch.Tensor

    @property
    def nnz(self) -> int:
        return self.qkeys.numel()


def make(cfg: Config, device="cpu", with_values: bool = True) -> Workload:
    keys = table_keys(cfg, device)
    offsets, qkeys = batch(cfg, device)
    n_elems = int(sum(cfg.vocab[s] * cfg.dims[s] for s in range(cfg.n_slots)))
    values = w0_values(cfg, n_elems, device) if with_values else None
    return Workload(cfg, keys, offsets, qkeys, values, grad_out(cfg, device))
