"""bench.py's recorded DRAM traffic (profiles/kda_traffic.json) on CPU: each kernel's figure is
reported only while the digest of that kernel's own sources matches the one recorded with it."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_every_recorded_kernel_has_its_source_list():
    with open(os.path.join(ROOT, "profiles", "kda_traffic.json")) as f:
        rec = json.load(f)
    assert set(rec["kernels"]) <= set(bench.KERNEL_SOURCES)
    for name, entry in rec["kernels"].items():
        assert entry["dram_bytes_per_launch"] > 0 and len(entry["source_sha256"]) == 64, name
        for src in bench.KERNEL_SOURCES[name]:
            assert os.path.exists(os.path.join(ROOT, "gated_delta_rule_08_gb300", "csrc", src)), src


def test_a_changed_source_drops_only_its_own_kernels(monkeypatch):
    real = bench.source_digest
    fresh = bench.measured_traffic()
    # pretend kda_decode.cu changed: only the decode kernel's traffic may disappear
    monkeypatch.setattr(bench, "source_digest",
                        lambda names: "0" * 64 if "kda_decode.cu" in names else real(names))
    after = bench.measured_traffic()
    assert "kda_decode" not in after
    assert {k: v for k, v in fresh.items() if k != "kda_decode"} == after


def test_digest_depends_on_names_and_contents():
    a = bench.source_digest(("kda_decode.cu", "kda_device.cuh"))
    b = bench.source_digest(("kda_device.cuh", "kda_decode.cu"))
    c = bench.source_digest(("kda_decode.cu",))
    assert len({a, b, c}) == 3
