"""Host logic of bench.py that needs no GPU: reading the committed ncu summary
of the scoring kernel for the roofline's traffic figure."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SCORE_SRC = os.path.join(ROOT, "sparse_attention_indexer_launch_gb300", "csrc", "score.cu")


def _summary_fields():
    fields = {}
    for line in open(os.path.join(ROOT, "profiles", "score_kernel_cfg3.md")):
        if line.startswith("- ") and ": " in line:
            k, v = line[2:].split(": ", 1)
            fields[k.strip()] = v.strip().strip("`")
    return fields


def test_summary_has_the_fields_bench_reads():
    f = _summary_fields()
    assert "score.cu sha256[:16]" in f
    assert int(f["dram bytes per launch"].replace(",", "")) > 0


def test_traffic_follows_the_kernel_source(tmp_path):
    import hashlib
    f = _summary_fields()
    sha = hashlib.sha256(open(SCORE_SRC, "rb").read()).hexdigest()[:16]
    got = bench.profile_traffic(SCORE_SRC)
    if f["score.cu sha256[:16]"] == sha:
        assert got == int(f["dram bytes per launch"].replace(",", ""))
    else:
        assert got is None
    # any other source text: the counters no longer describe it
    other = tmp_path / "score.cu"
    other.write_bytes(open(SCORE_SRC, "rb").read() + b"\n// changed\n")
    assert bench.profile_traffic(str(other)) is None


def test_cpu_baseline_sample_is_bounded_and_described():
    import oracle
    import workloads
    prob = workloads.make_config(0)           # one row of 4,096 keys: the oracle takes milliseconds
    orc = oracle.default()
    r = bench.cpu_baseline(prob, orc, budget_s=0.3)
    assert r["kind"] == "oracle" and r["unit"] == "key·rows/s"
    assert r["value"] > 0 and r["cores"] >= 1
    assert r["seconds"] < 2.0                 # about the budget, never far past it
    assert "pass(es) over the whole workload" in r["sample"]   # the workload fits: whole passes
    # a budget far below one pass cuts the rows instead of repeating them
    cut = bench.cpu_baseline(prob, orc, budget_s=1e-7, rate_hint=r["rate"])
    assert "of 1 rows" in cut["sample"] and cut["value"] > 0
