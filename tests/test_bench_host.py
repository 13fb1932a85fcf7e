"""Host logic of bench.py that needs no GPU: the algorithmic byte and flop
counts behind the roofline, and the source-hash rule for recorded traffic."""
import hashlib
import json
import os

import pytest

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_resident_step_bytes(bench):
    """Every entry resident: the resolve reads and writes each 1152-byte row once
    (plus 12 bytes of ids per entry); the decode reads each row once, q, out, lse
    and 8 bytes of ids per entry; 151.8 MB and 84.95 MB per step."""
    w = W.WORKLOADS["resident"]
    n = w.B * w.K
    r_hbm, r_link, d_bytes, flops = bench.algorithmic(w, (n, 0, 0))
    assert r_hbm == n * 1152 * 2 + n * 12 and r_link == 0
    assert abs(r_hbm / 1e6 - 151.8) < 0.1
    q, out = w.B * w.H * 576 * 2, w.B * w.H * (512 * 2 + 4)
    assert d_bytes == n * 1152 + q + out + n * 8
    assert abs(d_bytes / 1e6 - 84.95) < 0.01
    assert flops == 2.0 * w.B * w.H * w.K * 1088


def test_misses_and_in_place(bench):
    w = W.WORKLOADS["noresident"]
    n, rb = w.B * w.K, w.row_bytes
    res, hot, miss = 0, n // 2, n - n // 2
    g = bench.algorithmic(w, (res, hot, miss))
    p = bench.algorithmic(w, (res, hot, miss), in_place=True)
    assert g[0] == hot * rb + n * rb + miss * rb + n * 12      # hits read, all written, slots
    assert p[0] == miss * rb + n * 12                          # only the slots
    assert g[1] == p[1] == miss * rb                            # host link: each miss once
    assert g[2] == p[2] and g[3] == p[3]                        # attention reads the same rows


def test_per_token_counts_distinct_rows_once(bench):
    """One list per query token: entries are B*T*K, but a row several tokens
    select is read once and a missing row crosses the link once."""
    w = W.WORKLOADS["hybrid"]
    entries = w.B * w.T * w.K
    distinct_rows, distinct_misses = 42606.0, 18320.0
    r_hbm, r_link, d_bytes, flops = bench.algorithmic(
        w, (500, 88000, 42000), in_place=True, per_token=(distinct_rows, distinct_misses))
    assert r_link == distinct_misses * w.row_bytes
    assert r_hbm == distinct_misses * w.row_bytes + entries * 12
    q, out = w.B * w.T * w.H * 576 * 2, w.B * w.T * w.H * (512 * 2 + 4)
    assert d_bytes == distinct_rows * w.row_bytes + q + out + entries * 8
    assert flops == 2.0 * w.B * w.T * w.H * w.K * 1088


def test_traffic_record_follows_the_source_hash(bench):
    """A recorded DRAM figure is reported only while the kernel's source is the
    one it was captured from, and only for the way rows reached attention in
    the capture (in place or gathered)."""
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for k in ("resolve", "decode"):
        src = rec[k]["source"]
        sha = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
        mode = rec[k]["in_place"]
        got = bench._traffic(k, src, mode)
        assert got == (rec[k]["dram_bytes_per_launch"] if sha == rec[k]["source_sha"] else None)
        assert bench._traffic(k, src, not mode) is None
