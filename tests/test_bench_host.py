"""Host-side logic of bench.py (CPU): the DRAM-traffic record of the roofline kernel."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def _record(tmp_path, sha, nbytes=1000, tokens=10):
    name, _ = bench.TRAFFIC_RECORDS["csa.attention"]
    (tmp_path / name).write_text(
        "# capture summary\n\n"
        f"- `traffic_bytes_per_launch`: `{nbytes}`\n"
        f"- `tokens_per_launch`: `{tokens}`\n"
        f"- `source_sha256`: `{sha}`\n")


def test_traffic_scaled_by_tokens_when_sources_match(tmp_path):
    sha = bench.kernel_source_hash(bench.TRAFFIC_RECORDS["csa.attention"][1])
    _record(tmp_path, sha, nbytes=1000, tokens=10)
    assert bench.measured_traffic("csa.attention", 80, str(tmp_path)) == 8000.0


def test_traffic_null_once_the_kernel_changed(tmp_path):
    _record(tmp_path, "0" * 64)
    assert bench.measured_traffic("csa.attention", 80, str(tmp_path)) is None


def test_traffic_null_without_a_record(tmp_path):
    assert bench.measured_traffic("csa.attention", 80, str(tmp_path)) is None
    assert bench.measured_traffic("hca.attention", 80) is None


def test_committed_record_parses():
    # the committed summary carries the three fields in the format the bench reads
    name, _ = bench.TRAFFIC_RECORDS["csa.attention"]
    text = open(os.path.join(os.path.dirname(bench.__file__), "profiles", name)).read()
    for key in ("traffic_bytes_per_launch", "tokens_per_launch", "source_sha256"):
        assert f"- `{key}`:" in text
