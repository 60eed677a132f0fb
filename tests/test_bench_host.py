"""Host-side logic of bench.py that needs no GPU: the lookup of captured DRAM traffic, which
the bench line may only report while the kernel's sources are the ones that were profiled."""
import hashlib
import json

import pytest

import bench


def _setup(root, src_text="kernel body v1\n", entries=None):
    (root / "profiles").mkdir()
    (root / "src").mkdir()
    src = root / "src" / "k.cu"
    src.write_text(src_text)
    digest = hashlib.sha256(src_text.encode()).hexdigest()
    if entries is None:
        entries = [{"kernel": "main_kernel", "workload": "w", "sources": {"src/k.cu": digest},
                    "dram_bytes_read": 1000, "dram_bytes_write": 24}]
    (root / "profiles" / "dram_traffic.json").write_text(json.dumps({"entries": entries}))
    return src


@pytest.fixture
def root(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_traffic_reported_while_sources_match(root):
    _setup(root)
    assert bench.captured_traffic("main_kernel", "w") == 1024


def test_traffic_stale_after_a_source_edit(root):
    src = _setup(root)
    src.write_text("kernel body v2\n")
    assert bench.captured_traffic("main_kernel", "w") is None


def test_traffic_stale_when_a_source_is_missing(root):
    src = _setup(root)
    src.unlink()
    assert bench.captured_traffic("main_kernel", "w") is None


def test_traffic_needs_the_same_kernel_and_workload(root):
    _setup(root)
    assert bench.captured_traffic("main_kernel", "other") is None
    assert bench.captured_traffic("other_kernel", "w") is None


def test_traffic_every_listed_source_must_match(root):
    src = _setup(root)
    second = root / "src" / "h.cuh"
    second.write_text("header\n")
    entries = [{"kernel": "main_kernel", "workload": "w",
                "sources": {"src/k.cu": hashlib.sha256(src.read_bytes()).hexdigest(),
                            "src/h.cuh": hashlib.sha256(b"older header\n").hexdigest()},
                "dram_bytes_read": 1, "dram_bytes_write": 1}]
    (root / "profiles" / "dram_traffic.json").write_text(json.dumps({"entries": entries}))
    assert bench.captured_traffic("main_kernel", "w") is None


def test_traffic_none_without_a_readable_file(root):
    assert bench.captured_traffic("main_kernel", "w") is None  # no profiles/ at all
    (root / "profiles").mkdir()
    (root / "profiles" / "dram_traffic.json").write_text("{ not json")
    assert bench.captured_traffic("main_kernel", "w") is None


def test_committed_entries_name_existing_sources_and_summaries():
    # every committed entry points at files of this repository and carries both byte counts
    import os
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        doc = json.load(f)
    assert doc["entries"]
    for e in doc["entries"]:
        assert e["dram_bytes_read"] > 0 and e["dram_bytes_write"] >= 0
        for rel in e["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, rel)), rel
        assert os.path.exists(os.path.join(bench.ROOT, e["summary"])), e["summary"]


def test_default_workload_dominant_kernel_traffic_is_current():
    # the default benchmark line reports the backward main kernel's DRAM traffic only while the
    # capture matches the committed sources: a kernel edit without a new capture fails here
    w = bench.W.WORKLOADS[5]
    kernel = "bwd_tc64_kernel" if w.d == 64 else "bwd_tc_kernel"
    assert bench.captured_traffic(kernel, w.name) is not None


def _clock_line(sm, mx=2070, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return f"0, {sm}, {mx}, 812.5, 0x0000000000000000, {hw}, {hwt}, {swt}, {cap}"


def test_clock_summary_median_and_no_reasons():
    c = bench.ClockSampler(0)
    c.lines = [_clock_line(2070), _clock_line(2055), _clock_line(2070)]
    c.first = 0
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}


def test_clock_summary_reports_throttle_reasons():
    c = bench.ClockSampler(0)
    c.lines = [_clock_line(1980, cap="Active"), _clock_line(1500, hwt="Active"), _clock_line(2070)]
    c.first = 0
    assert c.summary()["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_summary_counts_only_the_timed_region():
    # samples before the timed region are left out, except the last one before it began
    c = bench.ClockSampler(0)
    c.lines = [_clock_line(900, hw="Active"), _clock_line(1000), _clock_line(2070), _clock_line(2070)]
    c.first = 2
    s = c.summary()
    assert s["samples"] == 3 and s["reasons"] == [] and s["sm_mhz"] == 2070.0


def test_clock_summary_skips_unreadable_rows():
    c = bench.ClockSampler(0)
    c.lines = ["0, [N/A], [N/A], [N/A], 0x0, Not Active, Not Active, Not Active, Not Active", "garbage",
               _clock_line(2040)]
    c.first = 0
    s = c.summary()
    assert s["samples"] == 1 and s["sm_mhz"] == 2040.0
    empty = bench.ClockSampler(0)
    assert empty.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_oracle_sample_block_is_part_of_a_causal_workload():
    # the CPU baseline times the leading n x n block of long heads; for causal attention the
    # first n query rows see only the first n keys, so the block's O, LSE and dQ rows are the
    # workload's own
    import numpy as np
    from oracle import ref
    r = np.random.default_rng(5)
    N, n, d = 300, 128, 16
    q, k, v, do = (r.standard_normal((N, d)) for _ in range(4))
    O, L = ref.forward_head(q, k, v, 0.25, True, rows=np.arange(n))
    Ob, Lb = ref.forward_head(q[:n], k[:n], v[:n], 0.25, True)
    assert np.allclose(O, Ob, rtol=0, atol=1e-13) and np.allclose(L, Lb, rtol=0, atol=1e-13)
    dq = ref.backward_head(q, k, v, do, 0.25, True, q_rows=np.arange(n))[0]
    dqb = ref.backward_head(q[:n], k[:n], v[:n], do[:n], 0.25, True)[0]
    assert np.allclose(dq, dqb, rtol=0, atol=1e-12)


def test_oracle_sample_counts_the_block_flops():
    w = bench.W.WORKLOADS[5]
    el, fl, heads, n = bench.oracle_sample(w, 0.0, max_heads=1, inp=_tiny_inputs(w))
    assert n == bench.SAMPLE_ROWS and heads == 1
    assert fl == 4 * n * n * w.d * 3.5 / 2


def _tiny_inputs(w):
    # the sampler reads only the leading block of each head: a tensor that long is enough
    import torch
    n = bench.SAMPLE_ROWS
    return {x: torch.randn(1, 1, n, w.d, generator=torch.Generator().manual_seed(i)).to(torch.bfloat16)
            for i, x in enumerate(("q", "k", "v", "do"))}
