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


def test_reference_arm_runs_without_the_product_library():
    """The oracle arm builds its inputs on the host (the oracle's block-manager
    model and the seeded host generator): it never loads libpagedkv.so, and it
    needs no GPU."""
    import json
    import subprocess
    code = ("import sys, json; sys.argv = ['bench.py', '--impl', 'reference', '--workload', "
            "'tiny', '--steps', '1', '--warmup', '0']; sys.path.insert(0, %r); import bench; "
            "bench.main(); maps = open('/proc/self/maps').read(); "
            "print(json.dumps({'product': 'libpagedkv' in maps, "
            "'oracle': '_liboracle' in maps}))" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = r.stdout.strip().splitlines()
    line, libs = json.loads(lines[-2]), json.loads(lines[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert libs == {"product": False, "oracle": True}


def test_host_case_matches_the_block_manager_model_workload():
    """The oracle arm's tables hold every context token: ceil(ctx / B) blocks
    per sequence, all distinct within a sequence, and the shared-prefix
    workload's sequences of one group share their prompt's full blocks."""
    for name in ("tiny", "opt13b", "shared_prefix"):
        hc = bench.host_case(name)
        B = hc["B"]
        for s, t in enumerate(hc["tables"]):
            assert len(t) == -(-int(hc["ctx"][s]) // B) and len(set(t)) == len(t)
    hc = bench.host_case("shared_prefix")
    p_len, _ = bench.W.prompt_and_suffix_lens(hc["spec"])
    g = hc["spec"].extra["per_group"]
    for gi, p in enumerate(p_len):
        full = int(p) // hc["B"]
        heads = {tuple(hc["tables"][gi * g + c][:full]) for c in range(g)}
        assert len(heads) == 1
