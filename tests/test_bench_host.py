"""Host logic of bench.py that needs no GPU: the DRAM traffic figure of the
roofline object is taken from an ncu summary only while the kernel sources it
names still have the recorded sha256 prefixes."""
import hashlib
import os

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "paged_kv_cache_92_gb300", "csrc")


def _prefix(name, n=16):
    with open(os.path.join(CSRC, name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:n]


def test_traffic_is_read_while_the_sources_match(tmp_path):
    s = tmp_path / "summary.md"
    s.write_text("traffic_bytes_per_launch: 123456\n"
                 f"source_sha256_prefix: pa_device.cuh={_prefix('pa_device.cuh')} "
                 f"pa_decode_tc.cu={_prefix('pa_decode_tc.cu', 12)}\n")
    assert bench.profiled_traffic(str(s)) == 123456


def test_traffic_is_dropped_once_a_source_changed(tmp_path):
    stale = "0" * 16 if _prefix("pa_device.cuh") != "0" * 16 else "1" * 16
    s = tmp_path / "summary.md"
    s.write_text("traffic_bytes_per_launch: 123456\n"
                 f"source_sha256_prefix: pa_decode_tc.cu={_prefix('pa_decode_tc.cu')} "
                 f"pa_device.cuh={stale}\n")
    assert bench.profiled_traffic(str(s)) is None


def test_traffic_needs_both_records(tmp_path):
    s = tmp_path / "summary.md"
    s.write_text("traffic_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic(str(s)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md")) is None
