"""bench.py's host-side bookkeeping, without a GPU: the stored ncu traffic is
reported only for the CUDA sources it was measured on, and the kernel count
per step follows the sort's digit width."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import sparse_ctr_embedding_gb300 as E  # noqa: E402


def test_stored_traffic_requires_matching_sources(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    wl, per = next(iter(rec["workloads"].items()))
    kernel, value = next(iter(per.items()))
    monkeypatch.setattr(bench, "kernel_fingerprint", lambda: rec["fingerprint"])
    assert bench.stored_traffic(wl, kernel) == value
    assert bench.stored_traffic(wl, "no_such_kernel") is None
    monkeypatch.setattr(bench, "kernel_fingerprint", lambda: "0" * 64)
    assert bench.stored_traffic(wl, kernel) is None


def test_fingerprint_is_stable():
    fp = bench.kernel_fingerprint()
    assert len(fp) == 64 and fp == bench.kernel_fingerprint()


def test_fingerprint_ignores_comments_only():
    a = 'int f(int x) { return x + 1; }  // one\n/* two */\nconst char* s = "//not a comment";\n'
    b = '// header\nint f(int x) { return x + 1; }\n\nconst char* s = "//not a comment";  /* tail */\n'
    assert bench.strip_comments(a) == bench.strip_comments(b)
    assert "//not a comment" in bench.strip_comments(a)
    assert bench.strip_comments(a) != bench.strip_comments(a.replace("x + 1", "x + 2"))


def test_launches_per_step_follow_the_digit_width():
    # placement (6) + recording forward, 5 launches per radix pass, reduce, fixup, and from
    # 2^24 lookups the fold kernel; the backward sorts rows within a slot: the largest
    # slot's key count sets the passes
    big = 1 << 24
    assert bench.launches_per_step(1_562_500, E.EMB_SORT_DIGIT_BITS, nnz=big) == 7 + 3 * 5 + 3   # 21 bits, 3 passes
    assert bench.launches_per_step(1_562_500, E.EMB_SORT_DIGIT_BITS, nnz=big - 1) == 7 + 3 * 5 + 2
    assert bench.launches_per_step(16_383, E.EMB_SORT_DIGIT_BITS) == 7 + 2 * 5 + 2        # 14 bits, 2 passes
    assert bench.launches_per_step(16_384, E.EMB_SORT_DIGIT_BITS) == 7 + 3 * 5 + 2        # 15 bits, 3 passes
    assert bench.launches_per_step(100, 7) == 7 + 1 * 5 + 2
    # the dedupe forward: placement, expand, the sort, dedupe pooling; the backward skips its sort
    assert bench.launches_per_step(1_562_500, E.EMB_SORT_DIGIT_BITS, dedup=True, nnz=big) == 7 + 3 * 5 + 1 + 3
