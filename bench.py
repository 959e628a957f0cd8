#!/usr/bin/env python
"""Benchmark of the embedding step on GB300: forward (probe + gather + pool)
and backward (dedupe + segmented reduce + Adagrad) over one CSR batch of a
seeded synthetic workload, through the C ABI.

Default workload: the large configuration (64 slots, 100M keys, dim 128,
float16 weights + float32 accumulators, batch 131,072, Zipf(1.1) bag lengths
in [1, 256], Zipf(1.1) ids, 5% absent keys, mean pooling).  Its inputs are far
larger than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=5, help="workload 1..5")
    ap.add_argument("--wdtype", default=None, choices=["f32", "f16", "f16m"],
                    help="weight storage instead of the workload's own (f16m: f32 master rows + f16 copy)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--fwd", default="fused", choices=["fused", "dedup"],
                    help="forward: the fused lookup + pooling (default), or the within-batch dedupe forward "
                         "(pairs sorted first, each unique row read once; the backward then skips its sort)")
    ap.add_argument("--vocab-div", type=int, default=1, help="shrink keys per slot (profiling a small case)")
    ap.add_argument("--batch-div", type=int, default=1, help="shrink the batch (profiling a small case)")
    ap.add_argument("--cpu-samples", type=int, default=2048,
                    help="samples of the batch the CPU-baseline oracle runs (bounded sample)")
    ap.add_argument("--ref-samples", type=int, default=128, help="samples per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--pipeline-depth", type=int, default=2,
                    help="buffer sets of the e2e leg's batch pipeline (uploads run up to depth - 1 batches ahead)")
    return ap.parse_args()


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (string and character literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


# The sources of the step's kernels and of the table they read (the forward, the
# backward, the host table build and the shared device code): a stored ncu figure
# is tied to these.  The batch pipeline and the device table build are host-side
# orchestration the captured kernels do not depend on.
STEP_SOURCES = ("emb_bwd.cu", "emb_fwd.cu", "emb_internal.cuh", "emb_table.cu")


def kernel_fingerprint() -> str:
    """sha256 of the step kernels' sources and the C ABI header with comments removed: ties a
    stored ncu figure to the code it measured (an edit of comments alone keeps it)."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_ctr_embedding_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in STEP_SOURCES]
    for f in files + [os.path.join(ROOT, "include", "emb_gb300.h")]:
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()


def stored_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu capture (profiles/dram_traffic.json),
    or None when absent or taken on other kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("fingerprint") != kernel_fingerprint():
        return None
    return d.get("workloads", {}).get(workload, {}).get(kernel)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init(args):
    import torch
    import torch.distributed as dist

    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(ws, x: float) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def launches_per_step(max_slot_keys: int, digit_bits: int, dedup: bool = False, nnz: int = 0) -> int:
    """Kernels this library launches for one forward (recording, or with dedupe) + one recorded bwd call.
    The backward sorts rows within a slot, so the pass count follows the largest slot; the fold kernel
    runs from 2^24 lookups."""
    bits = max(1, int(max_slot_keys).bit_length())
    passes = max(1, math.ceil(bits / digit_bits))
    fold = 1 if nnz >= (1 << 24) else 0
    # placement (transpose + 3 scan kernels + region setup + tile map); recording fwd, or expand + the
    # sort + dedupe pooling; (count + 3 scan + scatter) per radix pass; reduce; fold; fixup
    if dedup:
        return 6 + 1 + passes * 5 + 1 + 2 + fold
    return 6 + 1 + passes * 5 + 2 + fold


# ------------------------------------------------------------------ oracle (CPU baseline / reference arm)

class OracleRunner:
    """The CPU oracle on bounded samples (prefixes of whole samples) of the batch."""

    def __init__(self, cfg, keys_np, off_np, q_np, grad_np):
        import numpy as np

        import oracle

        self.np = np
        self.oracle = oracle
        self.cfg = cfg
        t0 = time.time()
        self.T = oracle.Table(keys_np, cfg.capacity, cfg.dims)
        self.build_s = time.time() - t0
        self.keys = keys_np
        self.off, self.q, self.grad = off_np, q_np, grad_np
        self.eoff = self.T.elem_offsets() if not cfg.uniform_dim else None

    def prepare(self, b0: int, b1: int):
        """Inputs for samples [b0, b1): a CSR sub-batch and the initial rows it touches."""
        import torch

        import workload as W

        np, cfg = self.np, self.cfg
        S = cfg.n_slots
        o = self.off[b0 * S:b1 * S + 1]
        q = self.q[o[0]:o[-1]]
        off = o - o[0]
        grad = self.grad[b0:b1]
        _, rows = self.T.resolve(q)
        rows = np.unique(rows[rows >= 0])
        dims_rows = np.array(cfg.dims, dtype=np.int64)[self.keys[rows] >> 48]
        if cfg.uniform_dim:
            eoff = torch.arange(0, (self.keys.size + 1) * cfg.dims[0], cfg.dims[0], dtype=torch.int64)
        else:
            eoff = torch.from_numpy(self.eoff)
        vals = W.w0_rows(cfg, eoff, torch.from_numpy(rows), torch.from_numpy(dims_rows)).numpy()
        row_map = np.full(self.keys.size, -1, dtype=np.int64)
        starts = np.concatenate([[0], np.cumsum(dims_rows)[:-1]]).astype(np.int64)
        row_map[rows] = starts
        return off, q, grad, vals, row_map

    def step(self, prep):
        """One oracle step on the sample: forward, per-key gradients, Adagrad. Returns seconds."""
        np, cfg, oracle = self.np, self.cfg, self.oracle
        off, q, grad, vals, row_map = prep
        t0 = time.perf_counter()
        self.T.forward(off, q, cfg.pool, cfg.wdtype, vals, row_map=row_map)
        uk, rows, goff, G, _ = self.T.backward(off, q, cfg.pool, grad)
        idx = np.concatenate([np.arange(row_map[r], row_map[r] + (goff[i + 1] - goff[i]))
                              for i, r in enumerate(rows)]) if rows.size else np.zeros(0, np.int64)
        oracle.adagrad(G, vals[idx], np.full(idx.size, cfg.acc0, np.float32), cfg.lr, cfg.eps)
        return time.perf_counter() - t0


def host_arrays(wl):
    return (wl.keys.cpu().numpy(), wl.offsets.cpu().numpy(), wl.qkeys.cpu().numpy(), wl.grad.cpu().numpy())


def run_reference(args):
    """--impl reference: the CPU oracle, timed on the host cores, on samples of the same workload."""
    import torch

    import workload as W

    ws, rank, local = dist_init(args)
    if rank != 0:
        return
    cfg = W.config(args.config)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if dev == "cuda":
        torch.cuda.set_device(local)
    keys = W.table_keys(cfg, dev).cpu().numpy()
    off_t, q_t = W.batch(cfg, dev)
    grad = W.grad_out(cfg, dev).cpu().numpy()
    runner = OracleRunner(cfg, keys, off_t.cpu().numpy(), q_t.cpu().numpy(), grad)
    b = max(1, min(args.ref_samples, cfg.batch))
    times, lookups = [], []
    for k in range(args.warmup + args.steps):
        b0 = (k * b) % max(1, cfg.batch - b + 1)
        prep = runner.prepare(b0, b0 + b)
        t = runner.step(prep)
        if k >= args.warmup:
            times.append(t)
            lookups.append(prep[1].size)
    total_t = sum(times)
    v = sum(lookups) / total_t
    line = {"metric": "embedding lookups/s (fwd+bwd step)", "value": v, "unit": "lookups/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total_t / len(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "sample_samples_per_step": b},
            "cpu_baseline": {"value": v, "unit": "lookups/s", "cores": 1, "kind": "oracle",
                             "sample": f"{b} samples x {cfg.n_slots} slots per step, rotating through the batch; "
                                       f"single-threaded oracle, {os.cpu_count()} cores available; "
                                       f"table build {runner.build_s:.1f}s untimed"},
            "e2e": {"value": v, "unit": "lookups/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def run_ours(args):
    import numpy as np
    import torch

    import workload as W
    import sparse_ctr_embedding_gb300 as E

    ws, rank, local = dist_init(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    E.build() if rank == 0 else None
    barrier(ws)
    E.build()
    cfg = W.config(args.config)
    if args.vocab_div > 1 or args.batch_div > 1:
        cfg = W.scaled(cfg, args.vocab_div, args.batch_div)
    if args.wdtype and args.wdtype != cfg.wdtype:
        cfg = dataclasses.replace(cfg, wdtype=args.wdtype, name=f"{cfg.name}/{args.wdtype}")
    stream = torch.cuda.current_stream()

    # ---- workload (generated on the device, keys copied to the host for the table build)
    t0 = time.time()
    keys = W.table_keys(cfg, dev)
    offsets, qkeys = W.batch(cfg, dev)
    grad = W.grad_out(cfg, dev)
    n_elems = int(sum(cfg.vocab[s] * cfg.dims[s] for s in range(cfg.n_slots)))
    values = W.w0_values(cfg, n_elems, dev)
    keys_h = keys.cpu()
    torch.cuda.synchronize()
    t_gen = time.time() - t0
    # the table prepared on the GPU from device keys (layout identical to the
    # host preparation below; built once without weights to time the build)
    t0 = time.time()
    try:
        E.emb_table_create_device(cfg.dims, cfg.wdtype, keys, capacity=cfg.capacity, acc_init=cfg.acc0).close()
        t_create_dev = time.time() - t0
    except E.EmbError as e:
        t_create_dev = f"not built: {e.name}"
    torch.cuda.empty_cache()
    t0 = time.time()
    tbl = E.emb_table_create(cfg.dims, cfg.wdtype, keys_h, values=values, capacity=cfg.capacity,
                             acc_init=cfg.acc0)
    t_create = time.time() - t0
    del values, keys
    torch.cuda.empty_cache()
    st = tbl.stats
    nnz = qkeys.numel()
    n_bags = offsets.numel() - 1
    out = torch.empty((cfg.batch, cfg.sum_dims), dtype=torch.float32, device=dev)
    wsb = torch.empty(E.emb_bwd_workspace_size(tbl, n_bags, nnz), dtype=torch.uint8, device=dev)

    # ---- algorithmic bytes of one step (the bytes the method must move)
    wsz = 2 if cfg.wdtype in ("f16", "f16m") else 4   # bytes of a row element the forward gathers
    _, rows = E.emb_resolve(tbl, qkeys)
    hit = rows >= 0
    dims_t = torch.tensor(cfg.dims, dtype=torch.int64, device=dev)
    d_occ = dims_t[qkeys >> 48]
    n_hits = int(hit.sum())
    gather_bytes = int((d_occ * hit).sum()) * wsz
    del rows, hit, d_occ
    p_bar = st["sum_probe"] / max(1, st["n_keys"])
    io_bytes = 8 * nnz + 16 * nnz * p_bar + 4 * cfg.batch * cfg.sum_dims + 8 * (n_bags + 1)
    fwd_bytes = io_bytes + gather_bytes

    fwd = E.emb_lookup_fwd_dedup if args.fwd == "dedup" else E.emb_lookup_fwd_record
    fwd_name = ("forward with dedupe (expand + sort + dedup_pool_kernel)" if args.fwd == "dedup"
                else "fwd_pool_kernel")

    def step():
        # the forward records each occurrence's resolved row for the backward
        fwd(tbl, offsets, qkeys, cfg.pool, wsb, out=out)
        E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz, cfg.pool, grad, cfg.lr, cfg.eps, wsb)

    step()
    uk = torch.empty(nnz, dtype=torch.int64, device=dev)
    nu = torch.zeros(1, dtype=torch.int64, device=dev)
    E.emb_bwd_unique_keys(tbl, wsb, uk, nu)
    n_unique = int(nu.item())
    d_u = dims_t[uk[:n_unique] >> 48]
    # per updated element: weights and accumulator read and written; a master-copy
    # table updates the f32 master and writes the element's f16 copy
    rmw_bytes = int(d_u.sum()) * (2 * 4 + 8 + 2 if cfg.wdtype == "f16m" else 2 * wsz + 8)
    del uk, d_u
    # the backward's bytes: the cached 4-byte row id of every occurrence (what
    # replaces the re-read of its key and the re-probe), the offsets, grad_out,
    # and the read-modify-write of the hit rows
    bwd_bytes = 4 * nnz + 8 * (n_bags + 1) + 4 * cfg.batch * cfg.sum_dims + rmw_bytes
    # algorithmic bytes per launch of each kernel (sort and partial sums are overhead)
    kernel_bytes = {
        fwd_name: fwd_bytes,
        "segreduce_update_kernel": 4 * cfg.batch * cfg.sum_dims + rmw_bytes,
    }
    flags = E.emb_check_device_flag(tbl)

    for _ in range(max(0, args.warmup - 1)):
        step()
    torch.cuda.synchronize()
    barrier(ws)
    clocks = Clocks(local)
    clocks.start()
    K = args.steps
    # per step: start, forward done, the backward's phases, backward call done
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3 + len(E.BWD_PHASES))] for _ in range(K)]
    for e in ev:                      # torch creates the CUDA event on first record
        for x in e:
            x.record(stream)
    torch.cuda.synchronize()
    for k in range(K):
        ev[k][0].record(stream)
        fwd(tbl, offsets, qkeys, cfg.pool, wsb, out=out)
        ev[k][1].record(stream)
        E.emb_bwd_phase_events(tbl, ev[k][2:-1])
        E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz, cfg.pool, grad, cfg.lr, cfg.eps, wsb)
        ev[k][-1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    E.emb_bwd_phase_events(tbl, [])
    total_ms = ev[0][0].elapsed_time(ev[K - 1][-1])
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[-1]) for e in ev)
    phase_ms = {name: statistics.mean(e[1 + i].elapsed_time(e[2 + i]) for e in ev)
                for i, name in enumerate(E.BWD_PHASES)}
    total_ms = max_over_ranks(ws, total_ms)
    ms_step = total_ms / K
    flags |= E.emb_check_device_flag(tbl)
    kernel_ms = {fwd_name: fwd_ms,
                 "radix sort (count + scan + scatter kernels)": phase_ms["sort"],
                 "segreduce_update_kernel": phase_ms["reduce"], "fixup_kernel": phase_ms["fixup"]}

    # ---- end to end through the C ABI: every step's CSR batch and grad_out are
    # copied in from pinned host memory and its pooled output copied back.  The
    # copies run on two copy streams into double buffers, overlapped with the
    # neighbouring steps (a loader feeding batches), and the timed region runs
    # from the first upload to the last download.
    e2e = None
    if not args.no_e2e:
        off_h = offsets.cpu().pin_memory()
        q_h = qkeys.cpu().pin_memory()
        g_h = grad.cpu().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()  # downloads are serialised on one stream
        h2d = off_h.numel() * 8 + q_h.numel() * 8 + g_h.numel() * 4
        d2h = out_h.numel() * 4
        # the library's batch pipeline: uploads of the next batch (copy stream) and
        # the pooled output's download (second copy stream) overlap the step
        pipe = E.Pipeline(tbl, n_bags, nnz, depth=args.pipeline_depth, upload_grad=True, stream=stream)

        def run_e2e(n_steps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            tickets = [pipe.submit(off_h, q_h, g_h)]
            for i in range(n_steps):
                if i + 1 < n_steps:
                    tickets.append(pipe.submit(off_h, q_h, g_h))
                pipe.forward(tickets[i], cfg.pool, out_h=out_h)
                pipe.backward_adagrad(tickets[i], cfg.lr, cfg.eps)
            pipe.wait(tickets[-1])
            torch.cuda.synchronize()
            return (time.perf_counter() - t0) * 1e3

        run_e2e(2)
        barrier(ws)
        Ke = max(3, K)   # as many steps as the device-timed leg: fill and drain weigh less
        e2e_ms = max_over_ranks(ws, run_e2e(Ke)) / Ke
        pipe.close()
        e2e = {"value": ws * nnz / (e2e_ms * 1e-3), "unit": "lookups/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "pipeline_depth": args.pipeline_depth,
               "path": "emb_pipeline (C ABI): pinned host CSR batch + grad_out uploaded on the pipeline's copy "
                       "stream, recording forward + recorded backward on the compute stream, pooled output "
                       "downloaded on its second copy stream; host wall clock from the first upload to the "
                       "last download"}

    peak, peak_src = peaks()
    fwd_gbs = fwd_bytes / (fwd_ms * 1e-3) / 1e9
    bwd_gbs = bwd_bytes / (bwd_ms * 1e-3) / 1e9
    single = {k: v for k, v in kernel_ms.items() if k in kernel_bytes}
    dom = max(single, key=single.get)
    dom_gbs = kernel_bytes[dom] / (kernel_ms[dom] * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": dom, "achieved": dom_gbs, "peak": peak, "unit": "GB/s",
            "frac": dom_gbs / peak, "traffic": stored_traffic(cfg.name, dom), "peak_source": peak_src,
            "algorithmic_bytes_per_launch": kernel_bytes[dom], "ms_per_launch": kernel_ms[dom]}
    kernels = {k: {"ms": v, "share": v / ms_step,
                   **({"algorithmic_gbs": kernel_bytes[k] / (v * 1e-3) / 1e9,
                       "frac_of_peak": kernel_bytes[k] / (v * 1e-3) / 1e9 / peak} if k in kernel_bytes else {})}
               for k, v in kernel_ms.items()}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        keys_np, off_np, q_np, g_np = keys_h.numpy(), offsets.cpu().numpy(), qkeys.cpu().numpy(), grad.cpu().numpy()
        runner = OracleRunner(cfg, keys_np, off_np, q_np, g_np)
        b = max(1, min(args.cpu_samples, cfg.batch))
        prep = runner.prepare(0, b)
        t = runner.step(prep)
        cpu = {"value": prep[1].size / t, "unit": "lookups/s", "cores": 1, "kind": "oracle",
               "sample": f"first {b} of {cfg.batch} samples ({prep[1].size} lookups, all {cfg.n_slots} slots): "
                         f"forward + per-key gradients + Adagrad in {t:.1f}s on 1 of {os.cpu_count()} host cores; "
                         f"oracle table build {runner.build_s:.1f}s untimed"}

    line = {
        "metric": "embedding lookups/s (fwd+bwd step)", "value": ws * nnz / (ms_step * 1e-3), "unit": "lookups/s",
        "n_gpus": ws, "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": cfg.name, "keys": cfg.n_keys, "slots": cfg.n_slots, "dim": cfg.dims[0]
                   if cfg.uniform_dim else list(cfg.dims), "weights": cfg.wdtype, "batch": cfg.batch,
                   "bags": n_bags, "nnz": nnz, "hits": n_hits, "unique_keys": n_unique, "pool": cfg.pool,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas" if ws > 1 else "single"},
        "samples_per_s": ws * cfg.batch / (ms_step * 1e-3),
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_lookups_per_s": nnz / (fwd_ms * 1e-3),
        "fwd_algorithmic_gbs": fwd_gbs, "bwd_algorithmic_gbs": bwd_gbs,
        "fwd_frac_nominal_8tbs": fwd_gbs / NOMINAL_HBM_GBS, "bwd_frac_nominal_8tbs": bwd_gbs / NOMINAL_HBM_GBS,
        "roofline": roof,
        "kernels": kernels,
        "fwd_roofline": {"achieved": fwd_gbs, "frac": fwd_gbs / peak, "algorithmic_bytes": fwd_bytes},
        "bwd_roofline": {"achieved": bwd_gbs, "frac": bwd_gbs / peak, "algorithmic_bytes": bwd_bytes},
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": K * launches_per_step(st["max_slot_keys"], E.EMB_SORT_DIGIT_BITS, args.fwd == "dedup", nnz),
        "clocks": clk, "device_flags": flags,
        "setup_s": {"generate": t_gen, "table_create": t_create, "table_create_device": t_create_dev},
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    tbl.close()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
