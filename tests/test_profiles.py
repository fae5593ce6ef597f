"""The committed DRAM-traffic records the bench line reports (no GPU).

bench.py looks up the attention kernel's DRAM traffic per launch in
profiles/traffic.txt under a hash of the attention sources; an edit to those
sources that is not followed by a new capture leaves the bench line's
`traffic` null.  This keeps the records in step with the code.
"""
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_traffic_records_match_the_attention_sources():
    sha = bench.src_sha()
    for workload in ("bass_b8", "bass_b8_e4m3", "draft_bass_b8"):
        t = bench.traffic_record(sha, workload)
        assert t is not None, f"no traffic record for {workload} at attention source hash {sha}"
        assert 5e7 < t < 5e8, (workload, t)


def test_traffic_record_lines_are_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.txt")) as fh:
        for ln in fh:
            f = ln.split()
            assert len(f) == 4 and f[0] == "attention", ln
            assert len(f[2]) == 12 and int(f[2], 16) >= 0, ln
            assert int(f[3]) > 0, ln
