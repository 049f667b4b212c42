"""The benchmark's evidence records on CPU: a DRAM-traffic record counts only
while the kernels' sources still hash to the value it was captured on, and
every committed record is of a workload the benchmark knows, with a
plausible size."""
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from newton_schulz_06_gb300 import inputs as I  # noqa: E402


def test_committed_traffic_records_are_well_formed():
    recs = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    assert recs
    for key, ent in recs.items():
        kernel, workload = key.split("@")
        I.workload(workload)                       # a workload bench.py knows
        current = ent["source_sha"] == bench.source_sha(ent["source_files"])
        got = bench.traffic_for(kernel, workload)
        # reported exactly while current, never once a source has changed
        assert got == (ent["bytes_per_launch_full_workload"] if current else None), key
        assert 0 < ent["bytes_per_launch_full_workload"] < 2 * ent["algorithmic_bytes_per_launch"]


def test_traffic_record_goes_stale_when_a_source_changes(tmp_path, monkeypatch):
    # a copy of the repository's sources and records, with one kernel file
    # edited after the capture
    for d in ("profiles", os.path.join("newton_schulz_06_gb300", "csrc")):
        shutil.copytree(os.path.join(ROOT, d), tmp_path / d)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # as if just captured on these sources
    rec_path = tmp_path / "profiles" / "traffic.json"
    recs = json.loads(rec_path.read_text())
    ent = recs["ns2_kernel<3>@square_4096_bf16"]
    ent["source_sha"] = bench.source_sha(ent["source_files"])
    rec_path.write_text(json.dumps(recs))
    assert bench.traffic_for("ns2_kernel<3>", "square_4096_bf16") == \
        ent["bytes_per_launch_full_workload"]
    src = tmp_path / "newton_schulz_06_gb300" / "csrc" / "ns2_kernels.cu"
    src.write_text(src.read_text() + "\n// edited\n")
    assert bench.traffic_for("ns2_kernel<3>", "square_4096_bf16") is None
    assert bench.traffic_for("ns2_kernel<2>", "no_such_workload") is None
