"""bench.py's host-side reading of the committed ncu summaries (no GPU): a
roofline traffic figure is used only while the summary's kernel source digest
matches the sources, and a workload without a summary has none."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def committed_lines(name):
    kv = {}
    for line in open(os.path.join(ROOT, "profiles", name)):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            kv[k.strip()] = v.strip().strip("`")
    return kv


def test_traffic_follows_the_digest():
    for wl, prof, src in (("opt13b", None, None), ("short", None, None),
                          ("prefill", "paged_prefill_tc_prefill.md", bench.PREFILL_SOURCES)):
        kv = committed_lines(prof or "paged_decode_main_%s.md" % wl)
        digest = bench.kernel_source_digest(src) if src else bench.kernel_source_digest()
        t = bench.profiled_traffic(wl, prof, src)
        if kv["kernel_source_sha256_16"] == digest:
            assert t == float(kv["dram_bytes_per_launch_full_size"])
        else:
            assert t is None


def test_stale_digest_or_missing_summary_gives_none(monkeypatch):
    assert bench.profiled_traffic("tiny") is None
    monkeypatch.setattr(bench, "kernel_source_digest", lambda files=None: "0" * 16)
    assert bench.profiled_traffic("opt13b") is None
    assert bench.profiled_traffic("prefill", "paged_prefill_tc_prefill.md",
                                  bench.PREFILL_SOURCES) is None
